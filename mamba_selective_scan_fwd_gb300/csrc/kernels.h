// Kernel argument blocks and launchers (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "tma.cuh"

namespace ss {

struct FwdArgs {
    const void *u, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias;
    const float* h0;  // initial state [Bsz][Dch][N], or null (zero)
    void* y;
    float* last_state;
    int64_t Bsz, L, Dch, N;
    int softplus;
    int a_is_log;     // A holds A_log: the scan uses A = -exp(A_log)
    int dtype;        // 0 f32, 1 f16, 2 bf16
    // chunk summaries, per summary index (layout of FPlan): the end state from
    // a zero start [.][CH][N] and the chunk's sum of delta_eff [.][CH]
    float* ws_fsum;
    float* ws_fsd;
    // pre-gate readout y0 = sum_n h C + D u, f32 [Bsz][L][Dch], stored by the
    // saving and checkpoint passes for the backward's dz when z is given
    // (null: not stored)
    float* y0;
    // tiles staged by TMA through the kernel's tensor maps (else by per-thread
    // asynchronous copies), and the library's device status word, where a
    // kernel that gave up waiting for a copy leaves kDevWaitTimeout
    int use_tma;
    int* status;
};

// A[d, n] of the scan: the input itself, or -exp(A_log) in the A_log form.
__device__ __forceinline__ float scan_A(const FwdArgs& a, int64_t i) {
    const float v = a.A[i];
    return a.a_is_log ? -expf(v) : v;
}

struct BwdArgs {
    FwdArgs f;        // forward inputs; f.y / f.last_state unused
    const void* dy;
    const float* dlast;  // incoming gradient of last_state [Bsz][Dch][N], or null (zero)
    float *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *ddelta_bias;
    float* dh0;          // gradient of the initial state [Bsz][Dch][N], or null
    // reverse chunk summaries per summary index: the carry a chunk passes back
    // from a zero incoming adjoint [.][CH][N] and the chunk's sum of delta_eff [.][CH]
    float* ws_rsum;
    float* ws_rsd;
    const float* ws_ckpt;  // sub-chunk start states (layout of ckpt_bytes)
    const float* y0;       // the forward's pre-gate readout, f32 [Bsz][L][Dch]
    float* ws_bc;     // per-tile dB/dC partials: [2][tiles][Bsz][L][N]
    float* ws_dA;     // per-part dA partials: [q][CH][N]
    float* ws_dD;     // per-part dD partials: [q][CH]
    float* ws_db;     // per-part ddelta_bias partials: [q][CH]
};

// One decoding step in place on the state (ss_decode_step).
struct DecodeArgs {
    const void *u, *delta, *B, *C, *z;  // u, delta, z: io [Bsz, Dch]; B, C: io [Bsz, N]
    const float *A, *D, *delta_bias;
    float* state;                       // [Bsz][Dch][N], read and rewritten
    void* y;                            // io [Bsz, Dch]
    int64_t Bsz, Dch, N;
    int softplus, a_is_log, dtype;
};

// Workspace layout of the backward (byte offsets, each 256-aligned).
struct BwdLayout {
    size_t fsum, fsd, rsum, rsd, ckpt, bc, dA, dD, db, total;
};

constexpr int kModeY = 0, kModeSummary = 1, kModeCkpt = 2, kModeYSave = 3;

// Block layout shared by the forward and backward scans.  A lane holds S
// states of two adjacent channels (a channel pair), so every B / C value it
// reads from shared memory serves two channels.  For N >= 16 a block has two
// warps that split the states of every channel; within a warp G = NPW / S
// adjacent lanes share a channel pair, NPW = N / warps being the warp's
// states.  S is 4 where the warp holds at least four states (the backward
// keeps an 8-step window of the lane's 2 S states in registers: 64 floats),
// else all of them.  A block covers 2 * 32 / G channels (16 for N = 32, 32
// for N = 8 and 16, 64 for N <= 4) of one batch row and one time chunk.
__host__ __device__ constexpr int scan_warps(int64_t N) { return N >= 16 ? 2 : 1; }
__host__ __device__ constexpr int lane_states(int64_t N) {
    return N / scan_warps(N) >= 4 ? 4 : (int)(N / scan_warps(N));
}
__host__ __device__ constexpr int64_t channels_per_block(int64_t N) {
    return 2 * 32 / (N / scan_warps(N) / lane_states(N));
}

constexpr int kSub = 8;  // steps between saved states (the backward's recompute window)
constexpr int kFwdRows = 32;  // steps per forward tile

// Launch plan.  A unit is one (batch row, channel tile): unit u = b tiles_b +
// tile.  Units are grouped into at most two segments; a segment cuts the time
// axis of each of its units into K chunks of Lc steps (the last may be
// shorter), and every kernel launch covers one segment, one block per (unit,
// chunk).  Each (unit, chunk) is a part with an index q (segment order, then
// unit, then chunk) that places its parameter-gradient partials; the parts
// of chunked segments (K > 1) also have a summary index that places their
// chunk summaries.
struct Seg {
    int64_t u_lo, nu;  // units u_lo .. u_lo + nu
    int64_t K, Lc;     // chunks per unit and their length (a multiple of 32)
    int64_t q0;        // part of (u_lo, chunk 0); part (u, k) = q0 + (u - u_lo) K + k
    int64_t s0;        // summary index of (u_lo, chunk 0), likewise (K > 1 only)
};
struct FPlan {
    int64_t tiles_b;   // channel tiles (sizes the per-tile dB / dC partials)
    int64_t slots;     // saved-state slots per sequence: one per kSub steps of L rounded up to 32
    int nseg;
    Seg seg[2];
    int64_t parts;     // parts over all segments
    int64_t sparts;    // parts of the chunked segments (entries of the summary arrays)
    int64_t Kmax;      // the largest K
};

constexpr int64_t kSMs = 152;                  // SMs of a GB300
constexpr int64_t kTargetWarps = 8 * kSMs;     // 8 warps on every SM keep each one's pipes busy
constexpr int64_t kFwdMinChunk = 128;

// Bytes of chunk summaries (end state and sum of delta_eff per channel) that a
// split of a plan that needs none may add: within the 2 MiB scratch of the
// no-allocation forward, so that splitting never takes a problem out of it.
constexpr int64_t kSplitSummaryMax = 2 << 20;

// Forward declaration: blocks of one round (below).
inline int64_t round_blocks(int64_t N);

// Cost of cutting nunits units into K chunks of their L steps, in units of
// one round of full-length blocks: the rounds of chunk blocks, each 1 / K as
// long (a partial round counted whole), plus the chunk summaries, about 0.6 of
// a main pass for K - 1 of the K chunks.
inline double chunk_cost(int64_t nunits, int64_t K, int64_t rb) {
    return (double)ceil_div(nunits * K, rb) / (double)K +
           0.6 * (double)nunits / (double)rb * (double)(K - 1) / (double)K;
}

// Chunking of nunits units that fills the GPU: K time chunks when nunits
// blocks make less than one round, chosen by chunk_cost among the counts that
// fill at least one round (at most kcap; chunks of at least kFwdMinChunk
// steps; the cost is taken at the chunk length rounded up to 32 steps).
inline void chunking(int64_t nunits, int64_t L, int64_t N, int64_t& K, int64_t& Lc, int64_t kcap = 1ll << 40) {
    const int64_t rb = round_blocks(N);
    int64_t kmax = ceil_div(L, kFwdMinChunk);
    if (kmax > kcap) kmax = kcap;
    if (kmax < 1) kmax = 1;
    auto length = [&](int64_t k) {
        const int64_t lc = ceil_div(ceil_div(L, k), 32) * 32;
        return lc < 32 ? (int64_t)32 : lc;
    };
    K = 1;
    Lc = length(1);
    if (nunits <= 0 || nunits >= rb) return;
    const int64_t kmin = ceil_div(rb, nunits);
    double best = 0.0;
    bool have = false;
    for (int64_t k = kmin < kmax ? kmin : kmax; k <= kmax && k <= 3 * kmin; k++) {
        const int64_t lc = length(k), keff = ceil_div(L, lc);
        const double c = chunk_cost(nunits, keff, rb);
        if (!have || c < best - 1e-9) {
            best = c;
            have = true;
            K = keff;
            Lc = lc;
        }
    }
}

// Blocks of one round: kTargetWarps warps, 8 on every SM.  The scan kernels
// are built for 8 resident warps per SM (4 two-warp or 8 one-warp blocks:
// their register budget), so a round is also what one wave of the GPU holds.
inline int64_t round_blocks(int64_t N) { return kTargetWarps / scan_warps(N); }

// A pure function of the sizes (the same sizes always plan the same way).
// One segment chunked to fill the GPU; or, when the units already fill it, one
// block per unit -- except that a count of units that is not a whole number
// of rounds leaves a last partial round: its blocks run as a wave of their
// own on part of the GPU (each SM's throughput does not grow past 8 resident
// warps, and falls below it).  Those last units mod round units then form a
// second segment cut in time, so that every SM gets an equal share, when that
// costs less than the partial round (estimated as at least half a round; the
// chunk summaries of the second segment take about 0.6 of a main pass).
inline FPlan make_fplan(int64_t Bsz, int64_t L, int64_t Dch, int64_t N) {
    FPlan p;
    p.tiles_b = ceil_div(Dch, channels_per_block(N));
    p.slots = ceil_div(L, 32) * (32 / kSub);
    const int64_t units = Bsz * p.tiles_b;
    p.nseg = 1;
    p.seg[0].u_lo = 0;
    p.seg[0].nu = units;
    p.seg[0].q0 = 0;
    p.seg[0].s0 = 0;
    chunking(units, L, N, p.seg[0].K, p.seg[0].Lc);
    p.seg[1] = p.seg[0];
    const int64_t rb = round_blocks(N);
    const int64_t tail = units % rb, rounds = units / rb;
    if (p.seg[0].K == 1 && tail > 0 && rounds > 0) {
        int64_t Kt, Lct;
        const int64_t kcap = kSplitSummaryMax / (tail * channels_per_block(N) * (N + 1) * 4);
        chunking(tail, L, N, Kt, Lct, kcap);
        if (Kt > 1) {
            // costs in rounds: the tail's chunks (whole rounds of them) and its summaries
            const double split = chunk_cost(tail, Kt, rb);
            const double partial = (double)tail / (double)rb > 0.5 ? (double)tail / (double)rb : 0.5;
            if (split < partial) {
                p.nseg = 2;
                p.seg[0].nu = units - tail;
                p.seg[1].u_lo = units - tail;
                p.seg[1].nu = tail;
                p.seg[1].K = Kt;
                p.seg[1].Lc = Lct;
                p.seg[1].q0 = units - tail;
            }
        }
    }
    p.parts = 0;
    p.sparts = 0;
    p.Kmax = 1;
    for (int i = 0; i < p.nseg; i++) {
        p.seg[i].s0 = p.sparts;
        p.parts += p.seg[i].nu * p.seg[i].K;
        if (p.seg[i].K > 1) p.sparts += p.seg[i].nu * p.seg[i].K;
        if (p.seg[i].K > p.Kmax) p.Kmax = p.seg[i].K;
    }
    return p;
}

// Segment si of the plan, by value (selected field by field, so that a
// kernel parameter is never indexed at run time).
__host__ __device__ inline Seg seg_at(const FPlan& p, int si) {
    Seg s;
    s.u_lo = si ? p.seg[1].u_lo : p.seg[0].u_lo;
    s.nu = si ? p.seg[1].nu : p.seg[0].nu;
    s.K = si ? p.seg[1].K : p.seg[0].K;
    s.Lc = si ? p.seg[1].Lc : p.seg[0].Lc;
    s.q0 = si ? p.seg[1].q0 : p.seg[0].q0;
    s.s0 = si ? p.seg[1].s0 : p.seg[0].s0;
    return s;
}

// Segment holding unit u.
__host__ __device__ inline Seg seg_of(const FPlan& p, int64_t u) {
    return seg_at(p, (p.nseg > 1 && u >= p.seg[1].u_lo) ? 1 : 0);
}

// Whether any segment is cut into chunks (the chunk summaries are needed).
inline bool plan_chunked(const FPlan& p) { return p.Kmax > 1; }


// Measurement aid behind ss_profile_events: prof_mark records the next of
// the caller's events on `st` (nothing when none are set); every launcher
// marks before each kernel it launches, the entry point once after the last.
void prof_mark(cudaStream_t st);

// Launchers of one io type T (float, __half, __nv_bfloat16), defined in the
// per-io translation units.
template <typename T>
cudaError_t launch_fwd_io(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt,
                          const TmaMaps& maps);
template <typename T>
cudaError_t launch_bwd_io(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out, const TmaMaps& fmaps,
                          const TmaMaps& bmaps);

// ckpt: where the Y-mode forward also stores the states entering every kSub-th step (may be null).
// maps: the forward's tensor maps (boxes of kFwdRows steps), used when a.use_tma.
cudaError_t launch_fwd(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt, const TmaMaps& maps);
// ckpt_out: the checkpoint buffer to fill first, or null when a.ws_ckpt already
// holds the states saved by the forward.
// fmaps / bmaps: tensor maps of the forward (checkpoint pass) and of the backward
// (boxes of kSub steps), used when a.f.use_tma.
cudaError_t launch_bwd(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out, const TmaMaps& fmaps,
                       const TmaMaps& bmaps);

// Carry pass of time-cut segment si (K > 1) in the backward, between the reverse
// summaries and the main pass: it folds the summaries into the adjoint carry
// into the end of every chunk, in place over the summaries the main pass reads.
cudaError_t launch_bwd_carry(const BwdArgs& a, const FPlan& p, int si, cudaStream_t st);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

// Bytes of what the forward keeps for the backward (ss_fwd_save writes it
// into the caller's buffer; ss_bwd's checkpoint pass into its workspace):
// the state entering every kSub-th step of every (b, d) row, which the
// backward recomputes its windows from, then at ckpt_y0_offset the pre-gate
// readout y0 (f32 [Bsz][L][Dch]).  States layout: [b][channel tile][slot t /
// kSub][block of CH x N floats] (ckpt_block): the blocks of consecutive slots
// of a unit are contiguous, so that the backward copies two at a time.
// Within a block, lane l of warp w holds S states of its first channel at
// ckpt_slot(w, l, S, 0) and S of its second at ckpt_slot(w, l, S, 1) (the
// scan kernels' lane layout): the 32 lanes' runs of one channel of their pair
// are contiguous, so that a warp's 16-byte stores and loads of them are 512
// contiguous bytes (and free of shared-memory bank conflicts once staged).
inline size_t ckpt_y0_offset(const FPlan& p, int64_t Bsz, int64_t N) {
    return align_up((size_t)Bsz * p.tiles_b * channels_per_block(N) * p.slots * N * sizeof(float), 256);
}
inline size_t ckpt_bytes(const FPlan& p, int64_t Bsz, int64_t L, int64_t Dch, int64_t N) {
    return ckpt_y0_offset(p, Bsz, N) + (size_t)Bsz * L * Dch * sizeof(float);
}

// Float offset of the saved-state block of (batch row b, channel tile, slot).
__host__ __device__ inline int64_t ckpt_block(const FPlan& p, int64_t b, int64_t tile, int64_t slot, int64_t N) {
    return ((b * p.tiles_b + tile) * p.slots + slot) * (channels_per_block(N) * N);
}

// Float offset of lane's S saved states of channel e (0: the first of its
// pair, 1: the second) within a saved-state block.
__host__ __device__ constexpr int64_t ckpt_slot(int w, int lane, int S, int e) {
    return ((int64_t)(2 * w + e) * 32 + lane) * S;
}

// Bytes of the forward chunk summaries (0 when nothing is chunked): end
// states [sparts][CH][N], then the sums of delta_eff [sparts][CH] at the
// 256-aligned offset fsum_offset_sd.
inline size_t fsum_offset_sd(const FPlan& p, int64_t N) {
    return align_up((size_t)p.sparts * channels_per_block(N) * N * sizeof(float), 256);
}
inline size_t fsum_bytes(const FPlan& p, int64_t N) {
    if (!plan_chunked(p)) return 0;
    return fsum_offset_sd(p, N) + align_up((size_t)p.sparts * channels_per_block(N) * sizeof(float), 256);
}

// Workspace of the backward (byte offsets, each 256-aligned): forward and
// reverse chunk summaries (only when chunked), sub-chunk start states (unless
// the forward saved them), per channel-tile dB / dC partials, per-part
// dA / dD / ddelta_bias partials.
inline BwdLayout bwd_layout2(const FPlan& p, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, bool saved) {
    BwdLayout w;
    size_t off = 0;
    const size_t pc = (size_t)p.parts * channels_per_block(N);    // partials
    const size_t sc = (size_t)p.sparts * channels_per_block(N);   // summaries
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    const bool ch = plan_chunked(p);
    w.fsum = take(ch && !saved ? sc * N * sizeof(float) : 0);
    w.fsd = take(ch && !saved ? sc * sizeof(float) : 0);
    w.rsum = take(ch ? sc * N * sizeof(float) : 0);
    w.rsd = take(ch ? sc * sizeof(float) : 0);
    w.ckpt = take(saved ? 0 : ckpt_bytes(p, Bsz, L, Dch, N));
    w.bc = take(2 * (size_t)p.tiles_b * Bsz * L * N * sizeof(float));
    w.dA = take(pc * N * sizeof(float));
    w.dD = take(pc * sizeof(float));
    w.db = take(pc * sizeof(float));
    w.total = off;
    return w;
}

}  // namespace ss
