// Kernel argument blocks and launchers (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

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
    int dtype;        // 0 f32, 2 bf16
    float* ws_fsum;   // chunk summaries (P, H): [Bsz*Dch][K][N] float2
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
    float* ws_rsum;   // reverse chunk summaries (P, M): [Bsz*Dch][K][N] float2
    const float* ws_ckpt;  // sub-chunk start states, step-major: [K * Lc/kSub][Bsz*Dch][N]
    float* ws_bc;     // per-tile dB/dC partials: [2][tiles][Bsz][L][N]
    float* ws_dA;     // per-(b,k) dA partials: [Bsz][K][Dch][N]
    float* ws_dD;     // per-(b,k) dD partials: [Bsz][K][Dch]
    float* ws_db;     // per-(b,k) ddelta_bias partials: [Bsz][K][Dch]
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
    size_t fsum, rsum, ckpt, bc, dA, dD, db, total;
};

constexpr int kModeY = 0, kModeSummary = 1, kModeCkpt = 2, kModeYSave = 3;

// Block layout shared by the forward and backward scans.  A lane holds S
// states of two adjacent channels (a channel pair), so every B / C value it
// reads from shared memory serves two channels.  For N >= 16 a block has two
// warps that split the states of every channel; within a warp G = 2 adjacent
// lanes share a channel pair (one lane for N = 1).  A block therefore covers
// 2 * 32 / G channels (32, or 64 for N = 1) of one batch row and one time
// chunk.
__host__ __device__ constexpr int fwd_warps(int64_t N) { return N >= 16 ? 2 : 1; }
__host__ __device__ constexpr int64_t channels_per_block(int64_t N) { return N >= 2 ? 32 : 64; }

// Launch plan: one block per (batch, channel tile, time chunk).  The time
// chunking (K, Lc) is shared by every kernel of a call.
struct FPlan {
    int64_t tiles_b; // channel tiles (sizes the per-tile dB / dC partials)
    int64_t K;       // time chunks
    int64_t Lc;      // chunk length (multiple of 32); the last chunk may be shorter
};

constexpr int64_t kTargetWarps = 1216;  // 8 warps on each of 152 SMs
constexpr int64_t kFwdMinChunk = 128;

// A pure function of the sizes (the same sizes always chunk the same way).
inline FPlan make_fplan(int64_t Bsz, int64_t L, int64_t Dch, int64_t N) {
    FPlan p;
    p.tiles_b = ceil_div(Dch, channels_per_block(N));
    const int64_t warps = Bsz * p.tiles_b * fwd_warps(N);
    int64_t K = 1;
    if (warps > 0 && warps < kTargetWarps) K = ceil_div(kTargetWarps, warps);
    const int64_t kmax = ceil_div(L, kFwdMinChunk);
    if (K > kmax) K = kmax;
    if (K < 1) K = 1;
    p.Lc = ceil_div(ceil_div(L, K), 32) * 32;
    if (p.Lc < 32) p.Lc = 32;
    p.K = ceil_div(L, p.Lc);
    if (p.K < 1) p.K = 1;
    return p;
}

constexpr int kSub = 4;  // backward sub-chunk: steps whose states stay in registers (checkpoint interval)

// Measurement aid behind ss_profile_events: prof_mark records the next of
// the caller's events on `st` (nothing when none are set); every launcher
// marks before each kernel it launches, the entry point once after the last.
void prof_mark(cudaStream_t st);

// Launchers of one io type T (float, __half, __nv_bfloat16), defined in the
// per-io translation units.
template <typename T>
cudaError_t launch_fwd2_io(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt);
template <typename T>
cudaError_t launch_bwd2_io(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out);

// ckpt: where the Y-mode forward also stores the sub-chunk start states (may be null).
cudaError_t launch_fwd2(const FwdArgs& a, const FPlan& p, cudaStream_t st, int mode, float* ckpt);
// ckpt_out: the checkpoint buffer to fill first, or null when a.ws_ckpt already
// holds the states saved by the forward.
cudaError_t launch_bwd2(const BwdArgs& a, const FPlan& p, cudaStream_t st, float* ckpt_out);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

// Bytes of the sub-chunk start states of every (b, d) row: the checkpoints the
// backward recomputes from (ss_fwd_save writes them into the caller's buffer).
// Layout: [k (Lc / kSub) + j][b][channel tile][block of CH x N floats]; within
// a block, float ((w 2 + e) 32 + lane) S + s is state n0 + s of channel c0 + e
// of the lane (the scan kernels' lane layout), so that a warp's stores and
// loads of one channel parity are contiguous.
inline size_t ckpt_bytes(const FPlan& p, int64_t Bsz, int64_t Dch, int64_t N) {
    (void)Dch;
    return (size_t)Bsz * p.tiles_b * channels_per_block(N) * p.K * (p.Lc / kSub) * N * sizeof(float);
}

// Float offset of a lane's slot for channel parity e within a saved-state block.
__host__ __device__ constexpr int64_t ckpt_slot(int w, int e, int lane, int S) {
    return ((int64_t)(w * 2 + e) * 32 + lane) * S;
}

// Workspace of the backward (byte offsets, each 256-aligned): forward and
// reverse chunk summaries (only when chunked), sub-chunk start states (unless
// the forward saved them), per channel-tile dB / dC partials, per-(batch,
// chunk) dA / dD / ddelta_bias partials.
inline BwdLayout bwd_layout2(const FPlan& p, int64_t Bsz, int64_t L, int64_t Dch, int64_t N, bool saved) {
    BwdLayout w;
    size_t off = 0;
    const size_t rows = (size_t)(Bsz * Dch);
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    w.fsum = take(p.K > 1 && !saved ? rows * p.K * N * 2 * sizeof(float) : 0);
    w.rsum = take(p.K > 1 ? rows * p.K * N * 2 * sizeof(float) : 0);
    w.ckpt = take(saved ? 0 : ckpt_bytes(p, Bsz, Dch, N));
    w.bc = take(2 * (size_t)p.tiles_b * Bsz * L * N * sizeof(float));
    w.dA = take((size_t)Bsz * p.K * Dch * N * sizeof(float));
    w.dD = take((size_t)Bsz * p.K * Dch * sizeof(float));
    w.db = take((size_t)Bsz * p.K * Dch * sizeof(float));
    w.total = off;
    return w;
}

}  // namespace ss
