// Launch dispatch on the io type (the kernels of each io type live in their
// own translation unit: fwd_*.cu, bwd_*.cu), and the backward's kernels that
// do not depend on it: the carry pass of time-cut segments and the two
// reductions.
#include "common.cuh"
#include "kernels.h"
#include "simd.cuh"

namespace ss {

// mode kModeY: the forward (summaries of the chunked segments, then y and
// last_state), also storing the state entering every kSub-th step into ckpt
// and the pre-gate readout into a.y0 when ckpt is given; mode kModeCkpt:
// the same walk writing only those states and the pre-gate readout (used by
// the backward), no y.
cudaError_t launch_fwd(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt, const TmaMaps& maps) {
    if (a.dtype == 0) return launch_fwd_io<float>(a, p, st, mode, ckpt, maps);
    if (a.dtype == 1) return launch_fwd_io<__half>(a, p, st, mode, ckpt, maps);
    return launch_fwd_io<__nv_bfloat16>(a, p, st, mode, ckpt, maps);
}

__global__ void k_bwd_reduce_bc(BwdArgs a, FPlan p);
__global__ void k_bwd_reduce_params(BwdArgs a, FPlan p);

// The backward's scan kernels (io-typed), then the two reductions.
cudaError_t launch_bwd(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out, const TmaMaps& fmaps,
                       const TmaMaps& bmaps) {
    cudaError_t e;
    if (a.f.dtype == 0) e = launch_bwd_io<float>(a, p, st, ckpt_out, fmaps, bmaps);
    else if (a.f.dtype == 1) e = launch_bwd_io<__half>(a, p, st, ckpt_out, fmaps, bmaps);
    else e = launch_bwd_io<__nv_bfloat16>(a, p, st, ckpt_out, fmaps, bmaps);
    if (e != cudaSuccess) return e;
    const int64_t n_bc = 2 * a.f.Bsz * a.f.L * a.f.N / (a.f.N % 4 == 0 ? 4 : 1);  // threads
    prof_mark(st);
    k_bwd_reduce_bc<<<(unsigned)ceil_div(n_bc, 256), 256, 0, st>>>(a, p);
    const int64_t n_par = a.f.Dch * a.f.N;
    prof_mark(st);
    k_bwd_reduce_params<<<(unsigned)ceil_div(n_par, 256), 256, 0, st>>>(a, p);
    return cudaGetLastError();
}

// Carry pass of a time-cut segment in the backward (one thread per (unit,
// channel, state)): from the reverse chunk summaries it forms the adjoint
// carry into the end of every chunk, so that a main-pass block reads its
// carry instead of folding the summaries of all the unit's later chunks
// itself.  r_{K-1} = d(last_state) (zero without one) and r_{k-1} = P_k r_k +
// M_k for k = K-1 .. 1, with M_k the carry chunk k passes back from a zero
// incoming adjoint and P_k = exp2(A log2(e) * the chunk's sum of delta_eff):
// each step is the one the main pass would take, in the same order and
// arithmetic, so the results are the same bits.  r_{k-1}, the carry into the
// end of chunk k - 1, is written over M_k, which nothing reads after it.  The
// summaries of eight chunks are loaded before they are folded, so that a
// thread waits for memory once per eight chunks.
constexpr int kCarryBatch = 8;

__global__ void k_bwd_carry(BwdArgs a, FPlan p, int si) {
    const FwdArgs& f = a.f;
    const Seg sgm = seg_at(p, si);
    const int64_t N = f.N, CH = channels_per_block(N), Dch = f.Dch;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= sgm.nu * CH * N) return;
    const int64_t ul = e / (CH * N), c = (e / N) % CH, n = e % N;
    const int64_t unit = sgm.u_lo + ul, b = unit / p.tiles_b, d = (unit % p.tiles_b) * CH + c;
    const bool ok = d < Dch;  // channels past Dch: read as zero by the main pass
    const float A2 = ok ? scan_A(f, d * N + n) * kLog2eF : 0.f;
    float r = ok && a.dlast ? a.dlast[(b * Dch + d) * N + n] : 0.f;
    const int64_t s_first = sgm.s0 + ul * sgm.K;         // reverse summaries of chunks 1 .. K-1
    float* M = a.ws_rsum + (s_first * CH + c) * N + n;  // chunk j at M[j CH N]
    const float* sd = a.ws_rsd + s_first * CH + c;     // chunk j at sd[j CH]
    for (int64_t j0 = sgm.K - 1; j0 >= 1; j0 -= kCarryBatch) {
        float mv[kCarryBatch], sv[kCarryBatch];
#pragma unroll
        for (int i = 0; i < kCarryBatch; i++) {
            const int64_t j = j0 - i >= 1 ? j0 - i : 1;  // below chunk 1: read, not folded
            mv[i] = M[j * CH * N];
            sv[i] = sd[j * CH];
        }
#pragma unroll
        for (int i = 0; i < kCarryBatch; i++) {
            if (j0 - i >= 1) {
                r = fmaf(ex2a(A2 * sv[i]), r, mv[i]);
                M[(j0 - i) * CH * N] = r;  // the carry into the end of chunk j0 - i - 1
            }
        }
    }
}

cudaError_t launch_bwd_carry(const BwdArgs& a, const FPlan& p, int si, cudaStream_t st) {
    const int64_t n = p.seg[si].nu * channels_per_block(a.f.N) * a.f.N;
    prof_mark(st);
    k_bwd_carry<<<(unsigned)ceil_div(n, 256), 256, 0, st>>>(a, p, si);
    return cudaGetLastError();
}

// dB / dC: sum of the per-tile partials, tiles in ascending order.  A thread
// owns 4 consecutive outputs (16-byte streaming loads, 8 tiles in flight)
// when N is a multiple of 4, one output otherwise.
__global__ void k_bwd_reduce_bc(BwdArgs a, FPlan p) {
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

// dA / dD / ddelta_bias: sum over the parts of each channel -- batch rows
// ascending, and within a row the chunks of its unit ascending.  The parts are
// visited in batches of kPB whose loads are all issued before their sums (the
// order of the sums is unchanged), so a thread waits for memory once per
// batch rather than once per part.
__global__ void k_bwd_reduce_params(BwdArgs a, FPlan p) {
    const int64_t Dch = a.f.Dch, N = a.f.N, CH = channels_per_block(N), Bsz = a.f.Bsz;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= Dch * N) return;
    const int64_t d = e / N, n = e % N;
    const int64_t tile = d / CH, c = d % CH;
    constexpr int kPB = 8;
    float acc = 0.f, accD = 0.f, accb = 0.f;
    int64_t b = 0, k = 0;  // the next part: chunk k of batch row b's unit
    Seg sg = seg_of(p, tile);
    while (b < Bsz) {
        int64_t qv[kPB];
#pragma unroll
        for (int j = 0; j < kPB; j++) {
            qv[j] = -1;
            if (b < Bsz) {
                qv[j] = sg.q0 + (b * p.tiles_b + tile - sg.u_lo) * sg.K + k;
                if (++k == sg.K) {
                    k = 0;
                    if (++b < Bsz) sg = seg_of(p, b * p.tiles_b + tile);
                }
            }
        }
        float v[kPB], vD[kPB], vb[kPB];
#pragma unroll
        for (int j = 0; j < kPB; j++) {
            v[j] = vD[j] = vb[j] = 0.f;
            if (qv[j] >= 0) {
                v[j] = a.ws_dA[(qv[j] * CH + c) * N + n];
                if (n == 0) {
                    vD[j] = a.ws_dD[qv[j] * CH + c];
                    vb[j] = a.ws_db[qv[j] * CH + c];
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kPB; j++) {
            if (qv[j] >= 0) {
                acc += v[j];
                accD += vD[j];
                accb += vb[j];
            }
        }
    }
    // A_log form: dA_log = dA * A with A = -exp(A_log)
    a.dA[e] = a.f.a_is_log ? acc * scan_A(a.f, e) : acc;
    if (n == 0) {
        if (a.dD) a.dD[d] = accD;
        if (a.ddelta_bias) a.ddelta_bias[d] = accb;
    }
}

}  // namespace ss
