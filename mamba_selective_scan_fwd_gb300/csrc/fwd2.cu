// Forward selective scan (baracuda-kernels `selective_scan.rs`, module doc
// "Algorithm summary"):
//
//   delta_eff = softplus?(delta + bias);  a = exp(delta_eff * A[d,n]);
//   h = a * h + delta_eff * B[t,n] * u;   y = (sum_n h * C[t,n] + D * u) * silu(z)
//
// One block owns CH channels of one batch row and one time chunk.  For
// N >= 16 the block has two warps and they split the N states of every
// channel: warp w holds states [w N/2, (w+1) N/2), G = 2 adjacent lanes per
// channel, S = N/4 states per lane.  Twice the warps of one-warp blocks keep
// the scheduler fed while each warp waits on MUFU and shared-memory results.
// Work per 32-step tile:
//   prologue  thread (warp w, lane l) takes time step t0 + l for channels
//             [w CH/NW, (w+1) CH/NW): converts its part of the row of u,
//             delta, z (contiguous runs of the [B, L, D] tensors), computes
//             delta_eff, delta_eff * u, silu(z) and D * u once per (t, d) and
//             stages them in shared memory; warp 0 stages the B row of its
//             step, warp 1 the C row;
//   scan      lane = (channel, state group) walks the 32 steps with packed
//             f32x2 arithmetic (one MUFU ex2 per state per step) and writes
//             its partial readout per step;
//   epilogue  thread (w, l) sums the partial readouts of step t0 + l over
//             the lanes and warps of each of its channels, adds D * u,
//             applies the gate and stores its part of the row of y.
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

template <typename T, int N>
struct FCfg {
    static constexpr int NW = fwd_warps(N);         // warps per block (they split the states)
    static constexpr int NPW = N / NW;              // states per warp
    static constexpr int G = NPW >= 2 ? 2 : 1;      // lanes per channel
    static constexpr int S = NPW / G;               // states per lane
    static constexpr int CH = 32 / G;               // channels per block
    static constexpr int CPT = CH / NW;             // channels per prologue / epilogue thread
    static constexpr int ESZ = (int)sizeof(T);
    static constexpr int RW = CPT * ESZ / 4;        // 32-bit words of a thread's part of a tile row
    static constexpr int NB = N * ESZ;              // bytes of a B / C row
    static constexpr int NWd = NB >= 4 ? NB / 4 : 1;  // 32-bit words per B / C row
    static constexpr int NP = N + 4;                // padded shared row of B / C (floats)
    static constexpr int YP = G == 2 ? 34 : 33;     // padded shared row of partial readouts
    static_assert(CPT * ESZ >= 16 && (CPT * ESZ) % 16 == 0, "a thread's row part is whole 16-byte vectors");
    static_assert(CH == kChannelsPerBlock || N == 1, "channel tile of the plan");
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

// CNT consecutive elements of a [Bsz, L, Dch] io tensor at element offset
// off (channel c0): vector loads when the run is aligned and complete,
// element loads (zero-filled past Dch) otherwise.
template <typename T, int CNT, int RW>
__device__ __forceinline__ void load_run(const T* base, int64_t off, int64_t c0, int64_t Dch, bool fast,
                                         uint32_t (&w)[RW]) {
    if (fast) {
        load_words<CNT * (int)sizeof(T), RW>(base + off, w);
    } else {
#pragma unroll
        for (int i = 0; i < RW; i++) w[i] = 0u;
#pragma unroll
        for (int c = 0; c < CNT; c++) {
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

// Stage a B or C row (N io elements held as words) as N floats of a shared row.
template <typename T, int N, int NWd>
__device__ __forceinline__ void stage_row(float* dst, const uint32_t (&w)[NWd], bool valid) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int n = 0; n < N; n += 4)
            *reinterpret_cast<float4*>(dst + n) =
                valid ? make_float4(elem<T>(w, n), elem<T>(w, n + 1), elem<T>(w, n + 2), elem<T>(w, n + 3))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
#pragma unroll
        for (int n = 0; n < N; n++) dst[n] = valid ? elem<T>(w, n) : 0.f;
    }
}

template <typename T, int N, int MODE>
__global__ void __launch_bounds__(32 * fwd_warps(N)) k_fwd2(FwdArgs a, FPlan p, int64_t ntiles, int64_t k_lo,
                                                            int64_t k_hi, float* ckpt) {
    constexpr bool SUMMARY = MODE == kModeSummary;
    constexpr bool NOY = MODE == kModeSummary || MODE == kModeCkpt;  // no readout, gate or y
    constexpr bool SAVE = MODE == kModeYSave || MODE == kModeCkpt;   // store the sub-chunk start states
    using C = FCfg<T, N>;
    constexpr int NW = C::NW, NPW = C::NPW, S = C::S, G = C::G, CH = C::CH, CPT = C::CPT, RW = C::RW,
                  NWd = C::NWd, NP = C::NP, YP = C::YP;
    // per-(t, d) staging, rows padded by one element: conflict-free for the
    // row-parallel prologue / epilogue (thread = step) and the scan (lane = channel)
    __shared__ float2 sDU[kRow][CH + 1];  // (delta_eff, delta_eff * u)
    __shared__ float2 sGD[NOY ? 1 : kRow][CH + 1];  // (gate, D * u)
    __shared__ __align__(16) float sB[kRow][NP];
    __shared__ __align__(16) float sC[NOY ? 1 : kRow][NP];
    __shared__ __align__(16) float sY[NOY ? 1 : NW][NOY ? 1 : kRow][YP];  // partial readouts, lane fastest
    __shared__ float sBias[CH], sDv[CH];

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
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

    if (tid < CH) {
        const int64_t dc = d0 + tid < Dch ? d0 + tid : Dch - 1;
        sBias[tid] = a.delta_bias ? a.delta_bias[dc] : 0.f;
        sDv[tid] = a.D ? a.D[dc] : 0.f;
    }

    // scan-lane identity: channel ch, states n0 .. n0 + S of warp w
    const int ch = lane / G, g = lane % G;
    const bool ch_ok = d0 + ch < Dch;
    const int64_t d = ch_ok ? d0 + ch : Dch - 1;
    const int n0 = w * NPW + g * S;
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
    // saved states, step-major: [k * (Lc / kSub) + j][Bsz * Dch][N]
    const int64_t ck_stride = a.Bsz * Dch * N;
    float* ck_row = SAVE ? ckpt + (k * (p.Lc / kSub)) * ck_stride + row * N + n0 : nullptr;

    // prologue-thread identity: step t0 + lane, channels cp0 .. cp0 + CPT
    const int cp0 = w * CPT;
    // B / C rows: with two warps, warp 0 stages B and warp 1 C; one warp stages both
    constexpr bool LOADB_ALL = NW == 1;
    const bool loads_b = LOADB_ALL || w == 0;
    const bool loads_c = !NOY && (LOADB_ALL || w == 1);
    uint32_t ru[RW], rd[RW], rz[RW], rb[NWd], rc[LOADB_ALL ? NWd : 1];
    auto load_rows = [&](int64_t t) {
        if (t < t_end) {
            const int64_t off = (b * L + t) * Dch + d0 + cp0;
            load_run<T, CPT, RW>(delta, off, d0 + cp0, Dch, fast, rd);
            load_run<T, CPT, RW>(u, off, d0 + cp0, Dch, fast, ru);
            if (!NOY && z) load_run<T, CPT, RW>(z, off, d0 + cp0, Dch, fast, rz);
            if constexpr (LOADB_ALL) {
                load_words<C::NB, NWd>(Bm + (b * L + t) * N, rb);
                if (!NOY) load_words<C::NB, NWd>(Cm + (b * L + t) * N, rc);
            } else {
                if (loads_b || loads_c) load_words<C::NB, NWd>((loads_b ? Bm : Cm) + (b * L + t) * N, rb);
            }
        }
    };
    load_rows(t_begin + lane);
    __syncthreads();

    for (int64_t t0 = t_begin; t0 < t_end; t0 += kRow) {
        // ---- prologue: step t0 + lane, channels cp0 .. cp0 + CPT
        {
            const bool rv = t0 + lane < t_end;
#pragma unroll
            for (int c = 0; c < CPT; c++) {
                const int cc = cp0 + c;
                float dl = 0.f, dlu = 0.f;
                if (rv) {
                    const float x = elem<T>(rd, c) + sBias[cc];
                    dl = a.softplus ? softplus_fast(x) : x;
                    dlu = dl * elem<T>(ru, c);
                }
                sDU[lane][cc] = make_float2(dl, dlu);
                if (!NOY) {
                    float gate = 1.f;
                    if (z) {
                        const float zz = elem<T>(rz, c);
                        gate = zz * sigmoid_fast(zz);
                    }
                    sGD[lane][cc] = make_float2(gate, sDv[cc] * elem<T>(ru, c));
                }
            }
            if constexpr (LOADB_ALL) {
                stage_row<T, N, NWd>(&sB[lane][0], rb, rv);
                if (!NOY) stage_row<T, N, NWd>(&sC[lane][0], rc, rv);
            } else {
                if (loads_b) stage_row<T, N, NWd>(&sB[lane][0], rb, rv);
                else if (loads_c) stage_row<T, N, NWd>(&sC[lane][0], rb, rv);
            }
        }
        if (t0 + kRow < t_end) load_rows(t0 + kRow + lane);
        __syncthreads();

        // ---- scan: 32 steps of this lane's S states.  Steps past t_end (last
        // tile only) carry delta_eff = 0 and B = 0: the state stays unchanged.
        float* ck_t = SAVE ? ck_row + ((t0 - t_begin) / kSub) * ck_stride : nullptr;
#pragma unroll 8
        for (int i = 0; i < kRow; i++) {
            if (SAVE && (i % kSub) == 0) {
                float* dst = ck_t + (i / kSub) * ck_stride;
                if constexpr (S % 4 == 0) {
#pragma unroll
                    for (int s = 0; s < S; s += 4)
                        if (ch_ok) *reinterpret_cast<float4*>(dst + s) = make_float4(h[s], h[s + 1], h[s + 2], h[s + 3]);
                } else {
#pragma unroll
                    for (int s = 0; s < S; s++)
                        if (ch_ok) dst[s] = h[s];
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
                if (!NOY) sY[w][i][lane] = yacc.x + yacc.y;
            } else {
                const float da = ex2a(du.x * A2[0]);
                h[0] = fmaf(da, h[0], du.y * Bv[0]);
                if (SUMMARY) P[0] *= da;
                else if (!NOY) sY[w][i][lane] = Cv[0] * h[0];
            }
        }
        __syncthreads();

        // ---- epilogue: step t0 + lane, channels cp0 .. cp0 + CPT
        if (!NOY) {
            const int64_t t = t0 + lane;
            if (t < t_end) {
                float yv[CPT];
#pragma unroll
                for (int c = 0; c < CPT; c++) {
                    const int cc = cp0 + c;
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < NW; q++) {
                        if constexpr (G == 2) {
                            const float2 v = *reinterpret_cast<const float2*>(&sY[q][lane][cc * 2]);
                            acc += v.x + v.y;
                        } else {
                            acc += sY[q][lane][cc];
                        }
                    }
                    const float2 gd = sGD[lane][cc];
                    yv[c] = (acc + gd.y) * gd.x;
                }
                T* yrow = static_cast<T*>(a.y) + (b * L + t) * Dch + d0 + cp0;
                if (fast) {
                    uint32_t wv[RW];
                    if constexpr (sizeof(T) == 4) {
#pragma unroll
                        for (int c = 0; c < CPT; c++) wv[c] = __float_as_uint(yv[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < CPT; c += 2) wv[c >> 1] = pack_bf16x2(yv[c], yv[c + 1]);
                    }
#pragma unroll
                    for (int v = 0; v < RW / 4; v++)
                        reinterpret_cast<uint4*>(yrow)[v] =
                            make_uint4(wv[4 * v], wv[4 * v + 1], wv[4 * v + 2], wv[4 * v + 3]);
                } else {
#pragma unroll
                    for (int c = 0; c < CPT; c++)
                        if (d0 + cp0 + c < Dch) st(yrow + c, yv[c]);
                }
            }
        }
    }

    if (SAVE && ch_ok) {
        // sub-chunk slots past the last tile (short last chunk only): the state
        // no longer changes there, so they hold the final state and the whole
        // buffer is written
        const int64_t nsub = p.Lc / kSub;
        const int64_t tiles_len = ((t_end - t_begin + kRow - 1) / kRow) * kRow;
        for (int64_t jj = tiles_len / kSub; jj < nsub; jj++) {
            float* dst = ck_row + jj * ck_stride;
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
    } else if (MODE != kModeCkpt && k == p.K - 1 && a.last_state && ch_ok) {
#pragma unroll
        for (int s = 0; s < S; s++) a.last_state[row * N + n0 + s] = h[s];
    }
}

template <typename T, int N>
int64_t fwd_tiles(int64_t Dch) {
    return ceil_div(Dch, FCfg<T, N>::CH);
}

template <typename T, int N, int MODE>
void launch_fwd_mode(const FwdArgs& a, const FPlan& p, cudaStream_t st, int64_t k_lo, int64_t k_hi, float* ckpt) {
    const int64_t nt = fwd_tiles<T, N>(a.Dch);
    prof_mark(st);
    k_fwd2<T, N, MODE><<<(unsigned)(nt * a.Bsz * (k_hi - k_lo)), 32 * FCfg<T, N>::NW, 0, st>>>(a, p, nt, k_lo,
                                                                                                 k_hi, ckpt);
}

template <typename T, int N>
cudaError_t launch_fwd2_t(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt) {
    if (p.K > 1) launch_fwd_mode<T, N, kModeSummary>(a, p, st, 0, p.K - 1, nullptr);
    if (mode == kModeCkpt) {
        launch_fwd_mode<T, N, kModeCkpt>(a, p, st, 0, p.K, ckpt);
    } else if (ckpt) {
        launch_fwd_mode<T, N, kModeYSave>(a, p, st, 0, p.K, ckpt);
    } else {
        launch_fwd_mode<T, N, kModeY>(a, p, st, 0, p.K, nullptr);
    }
    return cudaGetLastError();
}

// mode kModeY: the forward (summaries when K > 1, then y and last_state),
// also storing the state at every kSub-step sub-chunk start into ckpt when
// ckpt is given; mode kModeCkpt: the same walk writing only those states
// (used by the backward), no y.
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
