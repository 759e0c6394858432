// Kernel argument blocks and launchers (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace ss {

struct FwdArgs {
    const void *u, *delta, *B, *C, *z;
    const float *A, *D, *delta_bias;
    void* y;
    float* last_state;
    int64_t Bsz, L, Dch, N;
    int softplus;
    int dtype;        // 0 f32, 2 bf16
    float* ws_fsum;   // chunk summaries (P, H): [Bsz*Dch][K][N] float2
};

struct BwdArgs {
    FwdArgs f;        // forward inputs; f.y / f.last_state unused
    const void* dy;
    float *du, *ddelta, *dA, *dB, *dC, *dD, *dz, *ddelta_bias;
    float* ws_rsum;   // reverse chunk summaries M: [Bsz*Dch][K][N]
    float* ws_ckpt;   // sub-chunk start states: [Bsz*Dch*G][K][nsub][S]
    float* ws_bc;     // per-tile dB/dC partials: [2][tiles][Bsz][L][N]
    float* ws_dA;     // per-(b,k) dA partials: [Bsz][K][Dch][N]
    float* ws_dD;     // per-(b,k) dD partials: [Bsz][K][Dch]
    float* ws_db;     // per-(b,k) ddelta_bias partials: [Bsz][K][Dch]
};

// Workspace layout of the backward (byte offsets, each 256-aligned).
struct BwdLayout {
    size_t fsum, rsum, ckpt, bc, dA, dD, db, total;
};

inline BwdLayout bwd_layout(const Plan& p, int64_t Bsz, int64_t L, int64_t Dch, int64_t N) {
    BwdLayout w;
    size_t off = 0;
    const size_t rows = (size_t)(Bsz * Dch);
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    w.fsum = take(p.K > 1 ? rows * p.K * N * 2 * sizeof(float) : 0);
    w.rsum = take(p.K > 1 ? rows * p.K * N * sizeof(float) : 0);
    w.ckpt = take(rows * p.K * p.nsub * N * sizeof(float));
    w.bc = take(2 * (size_t)p.tiles * Bsz * L * N * sizeof(float));
    w.dA = take((size_t)Bsz * p.K * Dch * N * sizeof(float));
    w.dD = take((size_t)Bsz * p.K * Dch * sizeof(float));
    w.db = take((size_t)Bsz * p.K * Dch * sizeof(float));
    w.total = off;
    return w;
}

cudaError_t launch_fwd(const FwdArgs& a, const Plan& p, cudaStream_t st);
cudaError_t launch_fwd_summary(const FwdArgs& a, const Plan& p, cudaStream_t st);
cudaError_t launch_bwd(const BwdArgs& a, const Plan& p, cudaStream_t st);

}  // namespace ss
