// Forward selective scan (baracuda-kernels `selective_scan.rs`, module doc
// "Algorithm summary"):
//
//   delta_eff = softplus?(delta + bias);  a = exp(delta_eff * A[d,n]);
//   h = a * h + delta_eff * B[t,n] * u;   y = (sum_n h * C[t,n] + D * u) * silu(z)
//
// One warp owns CH = 32 / G channels of one batch row and one time chunk.
// Work per 32-step tile:
//   prologue  lane l takes time step t0 + l for all CH channels: converts the
//             row of u, delta, z (one contiguous CH-element run of the
//             [B, L, D] tensors) and the B / C rows, computes delta_eff,
//             delta_eff * u, silu(z) and D * u once per (t, d), and stages
//             them in shared memory;
//   scan      lane = (channel, state group): G lanes share a channel, each
//             holding S = N / G states in registers, and walk the 32 steps
//             with packed f32x2 arithmetic (one MUFU ex2 per state per step);
//   epilogue  lane l sums the G partial readouts of step t0 + l, adds D * u,
//             applies the gate and stores the row of y.
// The next tile's rows are loaded into registers while the current one is
// scanned.  The time axis is cut into K chunks only when batch x channels
// cannot fill the GPU; a chunk summary (P, H) = (product of a, end state
// from zero) then gives the carry-in state of the chunks after it.
#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"

namespace ss {

constexpr int kRow = 32;  // time steps per tile
static_assert(kRow % kSub == 0, "a tile holds whole checkpoint sub-chunks");

template <typename T, int N, int MODE>
struct FCfg {
    static constexpr int S = fwd_states_per_lane(N, MODE);  // states per lane
    static constexpr int G = N / S;                 // lanes per channel
    static constexpr int CH = 32 / G;               // channels per warp
    static constexpr int ESZ = (int)sizeof(T);
    static constexpr int ROWB = CH * ESZ;           // bytes of a tile row of a [B, L, D] tensor
    static constexpr int RW = ROWB / 4;             // 32-bit words per tile row
    static constexpr int NB = N * ESZ;              // bytes of a B / C row
    static constexpr int NW = NB >= 4 ? NB / 4 : 1; // 32-bit words per B / C row
    static constexpr int NP = N + 4;                // padded shared row of B / C (floats)
    static constexpr int YP = 32 + 4;               // padded shared row of partial readouts
};

// element j of a row held as 32-bit words
template <typename T>
__device__ __forceinline__ float elem(const uint32_t* w, int j) {
    if constexpr (sizeof(T) == 4) {
        return __uint_as_float(w[j]);
    } else {
        return (j & 1) ? bf16hi(w[j >> 1]) : bf16lo(w[j >> 1]);
    }
}

// Load NBYTES contiguous bytes (naturally aligned) into words.
template <int NBYTES, int NWORDS>
__device__ __forceinline__ void load_words(const void* p, uint32_t (&w)[NWORDS]) {
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

// Tile row of a [Bsz, L, Dch] io tensor at (b, t, d0..d0+CH): vector loads
// when the row is aligned and complete, element loads (zero-filled past Dch)
// otherwise.
template <typename T, int CH, int RW>
__device__ __forceinline__ void load_tile_row(const T* base, int64_t off, int64_t d0, int64_t Dch, bool fast,
                                              uint32_t (&w)[RW]) {
    if (fast) {
        load_words<CH * (int)sizeof(T), RW>(base + off, w);
    } else {
#pragma unroll
        for (int i = 0; i < RW; i++) w[i] = 0u;
#pragma unroll
        for (int c = 0; c < CH; c++) {
            if (d0 + c < Dch) {
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

// S consecutive floats of a shared row; the start is a multiple of S floats
// from a 16-byte aligned row, so S = 4, 8 use 16-byte loads.
template <int S>
__device__ __forceinline__ void ld_shared_row(const float* p, float (&v)[S]) {
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

template <typename T, int N, int MODE>
__global__ void __launch_bounds__(32) k_fwd2(FwdArgs a, FPlan p, int64_t ntiles, int64_t k_lo, int64_t k_hi,
                                             float* ckpt) {
    constexpr bool SUMMARY = MODE == kModeSummary;
    constexpr bool CKPT = MODE == kModeCkpt;
    constexpr bool NOY = SUMMARY || CKPT;  // no readout, gate or y
    using C = FCfg<T, N, MODE>;
    constexpr int S = C::S, G = C::G, CH = C::CH, RW = C::RW, NW = C::NW, NP = C::NP, YP = C::YP;
    // per-(t, d) staging, rows padded by one element: conflict-free for the
    // row-parallel prologue / epilogue (lane = step) and the scan (lane = channel)
    __shared__ float2 sDU[kRow][CH + 1];  // (delta_eff, delta_eff * u)
    __shared__ float2 sGD[kRow][CH + 1];  // (gate, D * u)
    __shared__ __align__(16) float sB[kRow][NP];
    __shared__ __align__(16) float sC[kRow][NP];
    __shared__ __align__(16) float sY[kRow][YP];
    __shared__ float sBias[CH], sDv[CH];

    const int lane = threadIdx.x;
    int64_t blk = blockIdx.x;
    const int64_t tile = blk % ntiles;
    blk /= ntiles;
    const int64_t nk = k_hi - k_lo;
    const int64_t k = k_lo + blk % nk;
    const int64_t b = blk / nk;
    const int64_t L = a.L, Dch = a.Dch;
    const int64_t d0 = tile * CH;
    const bool fast = ((Dch * (int64_t)sizeof(T)) % 16 == 0) && (d0 + CH <= Dch);
    const T* u = static_cast<const T*>(a.u);
    const T* delta = static_cast<const T*>(a.delta);
    const T* Bm = static_cast<const T*>(a.B);
    const T* Cm = static_cast<const T*>(a.C);
    const T* z = static_cast<const T*>(a.z);

    if (lane < CH) {
        const int64_t dc = d0 + lane < Dch ? d0 + lane : Dch - 1;
        sBias[lane] = a.delta_bias ? a.delta_bias[dc] : 0.f;
        sDv[lane] = a.D ? a.D[dc] : 0.f;
    }

    // scan-lane identity
    const int ch = lane / G, g = lane % G;
    const bool ch_ok = d0 + ch < Dch;
    const int64_t d = ch_ok ? d0 + ch : Dch - 1;
    const int n0 = g * S;
    float A2[S], h[S], P[S];
#pragma unroll
    for (int s = 0; s < S; s++) {
        A2[s] = a.A[d * N + n0 + s] * kLog2eF;
        h[s] = 0.f;
        P[s] = 1.f;
    }
    const int64_t row = b * Dch + d;
    if (!SUMMARY && k > 0) {
        const float2* sm = reinterpret_cast<const float2*>(a.ws_fsum) + row * p.K * N + n0;
        for (int64_t j = 0; j < k; j++) {
#pragma unroll
            for (int s = 0; s < S; s++) {
                const float2 ph = sm[j * N + s];
                h[s] = fmaf(ph.x, h[s], ph.y);
            }
        }
    }

    const int64_t t_begin = k * p.Lc;
    const int64_t t_end = t_begin + p.Lc < L ? t_begin + p.Lc : L;

    uint32_t ru[RW], rd[RW], rz[RW], rb[NW], rc[NW];
    auto load_rows = [&](int64_t t) {
        if (t < t_end) {
            const int64_t off = (b * L + t) * Dch + d0;
            load_tile_row<T, CH, RW>(delta, off, d0, Dch, fast, rd);
            load_tile_row<T, CH, RW>(u, off, d0, Dch, fast, ru);
            if (!NOY && z) load_tile_row<T, CH, RW>(z, off, d0, Dch, fast, rz);
            load_words<C::NB, NW>(Bm + (b * L + t) * N, rb);
            if (!NOY) load_words<C::NB, NW>(Cm + (b * L + t) * N, rc);
        }
    };
    load_rows(t_begin + lane);
    __syncwarp();

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kRow) {
        // ---- prologue: step t0 + lane, all CH channels
        {
            const bool rv = t0 + lane < t_end;
#pragma unroll
            for (int c = 0; c < CH; c++) {
                float dl = 0.f, dlu = 0.f;
                if (rv) {
                    const float x = elem<T>(rd, c) + sBias[c];
                    dl = a.softplus ? softplus_fast(x) : x;
                    dlu = dl * elem<T>(ru, c);
                }
                sDU[lane][c] = make_float2(dl, dlu);
                if (!NOY) {
                    float gate = 1.f;
                    if (z) {
                        const float zz = elem<T>(rz, c);
                        gate = zz * sigmoid_fast(zz);
                    }
                    sGD[lane][c] = make_float2(gate, sDv[c] * elem<T>(ru, c));
                }
            }
#pragma unroll
            for (int n = 0; n < N; n++) {
                sB[lane][n] = rv ? elem<T>(rb, n) : 0.f;
                if (!NOY) sC[lane][n] = rv ? elem<T>(rc, n) : 0.f;
            }
        }
        if (t0 + kRow < t_end) load_rows(t0 + kRow + lane);
        __syncwarp();

        // ---- scan: 32 steps of this lane's S states
#pragma unroll 8
        for (int i = 0; i < kRow; i++) {
            if (ckpt && (i % kSub) == 0 && ch_ok && t0 + i < t_end) {
                // state at the start of sub-chunk j = (t0 + i - t_begin) / kSub of chunk k,
                // stored step-major: [k * (Lc / kSub) + j][Bsz * Dch][N]
                const int64_t j = k * (p.Lc / kSub) + (t0 + i - t_begin) / kSub;
                float* dst = ckpt + (j * a.Bsz * a.Dch + row) * N + n0;
                if constexpr (S % 4 == 0) {
#pragma unroll
                    for (int s = 0; s < S; s += 4)
                        *reinterpret_cast<float4*>(dst + s) = make_float4(h[s], h[s + 1], h[s + 2], h[s + 3]);
                } else {
#pragma unroll
                    for (int s = 0; s < S; s++) dst[s] = h[s];
                }
            }
            const float2 du = sDU[i][ch];
            float Bv[S], Cv[S];
            ld_shared_row<S>(&sB[i][n0], Bv);
            if (!NOY) ld_shared_row<S>(&sC[i][n0], Cv);
            if constexpr (S >= 2) {
                const float2 dl2 = splat2(du.x), dlu2 = splat2(du.y);
                float2 yacc = make_float2(0.f, 0.f);
#pragma unroll
                for (int s = 0; s < S; s += 2) {
                    const float2 e = mul2(dl2, make_float2(A2[s], A2[s + 1]));
                    const float2 da = make_float2(ex2a(e.x), ex2a(e.y));
                    const float2 x = mul2(dlu2, make_float2(Bv[s], Bv[s + 1]));
                    const float2 hh = fma2(da, make_float2(h[s], h[s + 1]), x);
                    h[s] = hh.x;
                    h[s + 1] = hh.y;
                    if (SUMMARY) {
                        const float2 pp = mul2(make_float2(P[s], P[s + 1]), da);
                        P[s] = pp.x;
                        P[s + 1] = pp.y;
                    } else if (!NOY) {
                        yacc = fma2(make_float2(Cv[s], Cv[s + 1]), hh, yacc);
                    }
                }
                if (!NOY) sY[i][lane] = yacc.x + yacc.y;
            } else {
                const float da = ex2a(du.x * A2[0]);
                h[0] = fmaf(da, h[0], du.y * Bv[0]);
                if (SUMMARY) P[0] *= da;
                else if (!NOY) sY[i][lane] = Cv[0] * h[0];
            }
        }
        __syncwarp();

        // ---- epilogue: step t0 + lane, all CH channels
        if (!NOY) {
            const int64_t t = t0 + lane;
            if (t < t_end) {
                float yv[CH];
#pragma unroll
                for (int c = 0; c < CH; c++) {
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < G; q++) acc += sY[lane][c * G + q];
                    const float2 gd = sGD[lane][c];
                    yv[c] = (acc + gd.y) * gd.x;
                }
                T* yrow = static_cast<T*>(a.y) + (b * L + t) * Dch + d0;
                if (fast) {
                    uint32_t w[RW];
                    if constexpr (sizeof(T) == 4) {
#pragma unroll
                        for (int c = 0; c < CH; c++) w[c] = __float_as_uint(yv[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < CH; c += 2) w[c >> 1] = pack_bf16x2(yv[c], yv[c + 1]);
                    }
#pragma unroll
                    for (int v = 0; v < RW / 4; v++)
                        reinterpret_cast<uint4*>(yrow)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < CH; c++)
                        if (d0 + c < Dch) st(yrow + c, yv[c]);
                }
            }
        }
    }

    if (ckpt && ch_ok) {
        // sub-chunk slots past the end of the sequence (short last chunk only):
        // the state no longer changes there, so they hold the final state and
        // the whole checkpoint buffer is written
        const int64_t nsub = p.Lc / kSub;
        for (int64_t jj = (t_end - t_begin + kSub - 1) / kSub; jj < nsub; jj++) {
            float* dst = ckpt + ((k * nsub + jj) * a.Bsz * a.Dch + row) * N + n0;
#pragma unroll
            for (int s = 0; s < S; s++) dst[s] = h[s];
        }
    }

    if (SUMMARY) {
        if (ch_ok) {
            float2* out = reinterpret_cast<float2*>(a.ws_fsum) + (row * p.K + k) * N + n0;
#pragma unroll
            for (int s = 0; s < S; s++) out[s] = make_float2(P[s], h[s]);
        }
    } else if (!CKPT && k == p.K - 1 && a.last_state && ch_ok) {
#pragma unroll
        for (int s = 0; s < S; s++) a.last_state[row * N + n0 + s] = h[s];
    }
}

template <typename T, int N, int MODE>
int64_t fwd_tiles(int64_t Dch) {
    return ceil_div(Dch, FCfg<T, N, MODE>::CH);
}

template <typename T, int N>
cudaError_t launch_fwd2_t(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt) {
    if (p.K > 1) {
        const int64_t nt = fwd_tiles<T, N, kModeSummary>(a.Dch);
        prof_mark(st);
        k_fwd2<T, N, kModeSummary><<<(unsigned)(nt * a.Bsz * (p.K - 1)), 32, 0, st>>>(a, p, nt, 0, p.K - 1, nullptr);
    }
    if (mode == kModeCkpt) {
        const int64_t nt = fwd_tiles<T, N, kModeCkpt>(a.Dch);
        prof_mark(st);
        k_fwd2<T, N, kModeCkpt><<<(unsigned)(nt * a.Bsz * p.K), 32, 0, st>>>(a, p, nt, 0, p.K, ckpt);
    } else {
        const int64_t nt = fwd_tiles<T, N, kModeY>(a.Dch);
        prof_mark(st);
        k_fwd2<T, N, kModeY><<<(unsigned)(nt * a.Bsz * p.K), 32, 0, st>>>(a, p, nt, 0, p.K, ckpt);
    }
    return cudaGetLastError();
}

// mode kModeY: the forward (summaries when K > 1, then y and last_state);
// mode kModeCkpt: the same walk writing the state at every kSub-step
// sub-chunk start into ckpt (used by the backward), no y.
cudaError_t launch_fwd2(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt) {
#define SS_FWD2_N(T)                                                  \
    switch (a.N) {                                                    \
        case 1: return launch_fwd2_t<T, 1>(a, p, st, mode, ckpt);     \
        case 2: return launch_fwd2_t<T, 2>(a, p, st, mode, ckpt);     \
        case 4: return launch_fwd2_t<T, 4>(a, p, st, mode, ckpt);     \
        case 8: return launch_fwd2_t<T, 8>(a, p, st, mode, ckpt);     \
        case 16: return launch_fwd2_t<T, 16>(a, p, st, mode, ckpt);   \
        case 32: return launch_fwd2_t<T, 32>(a, p, st, mode, ckpt);   \
        default: return cudaErrorInvalidValue;                        \
    }
    if (a.dtype == 0) { SS_FWD2_N(float) }
    SS_FWD2_N(__nv_bfloat16)
#undef SS_FWD2_N
}

}  // namespace ss
